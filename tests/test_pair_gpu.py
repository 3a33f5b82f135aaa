"""Parity of the CTA-pair prefill kernel (FA_FLAG_PAIR: two-CTA clusters,
256-row MMAs, each CTA loading half of every K/V tile) with the fp64 oracle,
through the C ABI.  Gate: oracle/gate.py."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_and_check, run_kernel, sample_rows

pytestmark = pytest.mark.gpu

PAIR = fa.FA_FLAG_PAIR


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _assert(r):
    assert r.passed, str(r)


CASES = [  # B, H, Sq, Skv, dtype, causal
    (1, 1, 2, 2, "bf16", True),        # one pair item, almost all rows padding
    (1, 2, 129, 129, "bf16", True),    # ragged, stage 1 empty
    (1, 1, 257, 257, "fp16", False),   # stage 1 starts in the follower's half
    (1, 1, 513, 513, "bf16", True),    # two pair items, the second one row
    (2, 3, 1000, 1000, "bf16", True),
    (1, 1, 100, 300, "fp16", True),    # Sq < Skv (bottom-right diagonal)
    (1, 1, 300, 100, "bf16", True),    # Sq > Skv: rows without a visible key
    (1, 1, 600, 129, "fp16", True),
    (2, 8, 1024, 1024, "bf16", False),
    (2, 8, 1024, 1024, "bf16", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_pair_edge_shapes(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 128, dt, causal, 21, qk_mult=2.0, flags=PAIR))


# more pair items than pairs: every cluster takes several items in turn
PERSISTENT = [
    (4, 48, 600, 129, "bf16", True),
    (8, 32, 300, 300, "bf16", False),
    (1, 64, 1024, 128, "fp16", True),
]


@pytest.mark.parametrize("case", PERSISTENT, ids=lambda c: "x".join(map(str, c)))
def test_pair_persistent_item_sequences(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 128, dt, causal, 22, flags=PAIR))


def test_pair_headline_sampled_rows():
    w = inputs.HEADLINE
    rows = sample_rows(w.B, w.H, w.Sq, per_head=8, extra=256, seed=4)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=PAIR))


def test_pair_long_causal_sampled_rows():
    w = inputs.LONG16K
    rows = sample_rows(w.B, w.H, w.Sq, per_head=24, extra=128, seed=5)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=PAIR))


def test_pair_repeat_and_switches_bitwise_identical():
    q, k, v = inputs.make_qkv(2, 4, 1500, 1500, 128, "bf16", 23, 4.0)
    o1, l1 = run_kernel(q, k, v, True, flags=PAIR)
    o2, l2 = run_kernel(q, k, v, True, flags=PAIR)
    o3, l3 = run_kernel(q, k, v, True, flags=PAIR | fa.FA_FLAG_NO_LPT)
    o4, l4 = run_kernel(q, k, v, True, flags=PAIR | fa.FA_FLAG_ALWAYS_RESCALE)
    for o, l in ((o2, l2), (o3, l3), (o4, l4)):
        assert torch.equal(o, o1) and torch.equal(l, l1)


def test_single_cta_flag_on_a_pair_by_default_shape():
    """The headline shape runs on pairs by default; FA_FLAG_SINGLE_CTA runs
    the single-CTA kernel, which passes the same gate."""
    w = inputs.HEADLINE
    rows = sample_rows(w.B, w.H, w.Sq, per_head=4, extra=128, seed=6)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=fa.FA_FLAG_SINGLE_CTA))


def test_pair_flag_ignored_where_it_does_not_apply():
    """D=64 and an explicit key split run the single-CTA kernel."""
    _assert(run_and_check(1, 2, 300, 300, 64, "bf16", True, 24, flags=PAIR))
    q, k, v = inputs.make_qkv(1, 2, 256, 2048, 128, "bf16", 25)
    need = fa.fa_workspace_bytes(1, 2, 256, 2048, 128, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = run_kernel(q, k, v, True, flags=PAIR, num_splits=4, workspace=ws)
    _assert(check(q, k, v, o, lse, True, "bf16"))


def test_pair_watchdog_reports_timeout_and_context_survives():
    q, k, v = inputs.make_qkv(1, 2, 512, 512, 128, "bf16", 26)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)
    try:
        fa.fa_fwd_ex(dq, dk, dv, flags=PAIR | fa.FA_FLAG_TEST_STALL)
        assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_device_status() == fa.FA_OK
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = run_kernel(q, k, v, False, flags=PAIR)
    _assert(check(q, k, v, o, lse, False, "bf16"))


def test_pair_exact_running_max_mode():
    """FA_FLAG_EXACT_MAX on pairs passes the gate, and rescaling on every
    tile changes no bit."""
    w = inputs.C2_X4_CAUSAL
    q, k, v = w.make()
    o1, l1 = run_kernel(q, k, v, w.causal, flags=PAIR | fa.FA_FLAG_EXACT_MAX)
    _assert(check(q, k, v, o1, l1, w.causal, w.dtype))
    o2, l2 = run_kernel(q, k, v, w.causal,
                        flags=PAIR | fa.FA_FLAG_EXACT_MAX | fa.FA_FLAG_ALWAYS_RESCALE)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_pair_concurrent_streams_bitwise_identical():
    q, k, v = inputs.make_qkv(2, 8, 1024, 1024, 128, "bf16", 27)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ref, lref = fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=PAIR)
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for s in streams:
        with torch.cuda.stream(s):
            outs.append(fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=PAIR, stream=s))
    torch.cuda.synchronize()
    for o, l in outs:
        assert torch.equal(o, ref) and torch.equal(l, lref)
    assert fa.fa_get_device_status() == fa.FA_OK


def test_pair_scheduler_slots_wrap_around():
    """1100 pair launches (more than the 1024 scheduler slots), interleaved
    with single-CTA launches that share the slots: every launch claims every
    item."""
    q, k, v = inputs.make_qkv(2, 32, 1024, 512, 128, "bf16", 28)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ref, lref = fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=PAIR)
    o, lse = torch.empty_like(ref), torch.empty_like(lref)
    for i in range(1100):
        if i % 100 == 99:
            o.zero_()
            lse.fill_(float("nan"))
        fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=PAIR, out=o, lse=lse)
        if i % 7 == 3:
            fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=fa.FA_FLAG_SINGLE_CTA)
        if i % 100 == 99:
            torch.cuda.synchronize()
            assert torch.equal(o, ref) and torch.equal(lse, lref), i
    assert fa.fa_get_device_status() == fa.FA_OK


@pytest.mark.parametrize("case", [(4, 16, 4096, 4096, False), (2, 32, 2048, 2048, True),
                                  (8, 16, 1000, 1000, True)],
                         ids=lambda c: "x".join(map(str, c)))
def test_pair_many_items_per_cta_match_single_cta_bitwise(case):
    """Many items per pair (the item ring wraps dozens of times) give the
    same bits as the single-CTA kernel, which computes every element in the
    same order.  The pair kernel frees an item-ring slot with a relaxed
    cluster arrive, ordered after the read of the slot only by its control
    dependency on the value read; a slot overwritten before a taker read it
    would hand that taker another item and change the output here."""
    B, H, S, _, causal = case
    q, k, v = inputs.make_qkv(B, H, S, S, 128, "bf16", 71)
    ref = run_kernel(q, k, v, causal, flags=fa.FA_FLAG_SINGLE_CTA)
    for _ in range(3):
        o, lse = run_kernel(q, k, v, causal, flags=fa.FA_FLAG_PAIR)
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
