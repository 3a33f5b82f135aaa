"""Parity of the CTA-pair prefill kernel with 64-key score tiles and two
score buffers per stage (FA_FLAG_PAIR64) with the fp64 oracle, through the C
ABI.  Gate: oracle/gate.py."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_and_check, run_kernel, sample_rows

pytestmark = pytest.mark.gpu

P64 = fa.FA_FLAG_PAIR64


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _assert(r):
    assert r.passed, str(r)


CASES = [  # B, H, Sq, Skv, dtype, causal
    (1, 1, 2, 2, "bf16", True),        # one pair item, almost all rows padding
    (1, 1, 64, 64, "bf16", False),     # one key tile
    (1, 1, 65, 65, "fp16", True),      # a ragged second tile
    (1, 2, 129, 129, "bf16", True),    # stage 1 empty
    (1, 1, 257, 257, "fp16", False),   # stage 1 starts in the follower's half
    (1, 1, 513, 513, "bf16", True),    # two pair items, the second one row
    (2, 3, 1000, 1000, "bf16", True),
    (1, 1, 100, 300, "fp16", True),    # Sq < Skv (bottom-right diagonal)
    (1, 1, 300, 100, "bf16", True),    # Sq > Skv: rows without a visible key
    (1, 1, 600, 129, "fp16", True),
    (1, 1, 600, 40, "bf16", False),    # fewer keys than one tile
    (2, 8, 1024, 1024, "bf16", False),
    (2, 8, 1024, 1024, "bf16", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_pair64_edge_shapes(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 128, dt, causal, 31, qk_mult=2.0, flags=P64))


# more pair items than pairs: every cluster takes several items in turn
PERSISTENT = [
    (4, 48, 600, 129, "bf16", True),
    (8, 32, 300, 300, "bf16", False),
    (1, 64, 1024, 128, "fp16", True),
    (4, 16, 2048, 2048, "bf16", True),
]


@pytest.mark.parametrize("case", PERSISTENT, ids=lambda c: "x".join(map(str, c)))
def test_pair64_persistent_item_sequences(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 128, dt, causal, 32, flags=P64))


def test_pair64_headline_sampled_rows():
    w = inputs.HEADLINE
    rows = sample_rows(w.B, w.H, w.Sq, per_head=16, extra=256, seed=7)
    assert rows.size >= 512
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=P64))


def test_pair64_long_causal_sampled_rows():
    w = inputs.LONG32K
    rows = sample_rows(w.B, w.H, w.Sq, per_head=64, extra=256, seed=8)
    assert rows.size >= 512
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=P64))


def test_pair64_repeat_and_switches_bitwise_identical():
    """Repeats, the plain item order and rescaling on every tile give the
    same bits (many items per pair: the item ring wraps)."""
    q, k, v = inputs.make_qkv(4, 16, 1500, 1500, 128, "bf16", 33, 4.0)
    o1, l1 = run_kernel(q, k, v, True, flags=P64)
    o2, l2 = run_kernel(q, k, v, True, flags=P64)
    o3, l3 = run_kernel(q, k, v, True, flags=P64 | fa.FA_FLAG_NO_LPT)
    o4, l4 = run_kernel(q, k, v, True, flags=P64 | fa.FA_FLAG_ALWAYS_RESCALE)
    for o, l in ((o2, l2), (o3, l3), (o4, l4)):
        assert torch.equal(o, o1) and torch.equal(l, l1)


@pytest.mark.parametrize("scale", [1.0, 1e-3], ids=["sharp", "flat"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_pair64_extreme_scales(scale, causal):
    """A sharp softmax (the reference max moves, the rescale waits for the
    previous PV) and a nearly flat one; V scaled by 1/4 as in the other
    kernels' tests."""
    q, k, v = inputs.make_qkv(1, 4, 1500, 1500, 128, "bf16", 34)
    v = v * 0.25
    o, lse = run_kernel(q, k, v, causal, flags=P64, scale=scale)
    _assert(check(q, k, v, o, lse, causal, "bf16", scale=scale))


@pytest.mark.parametrize("exact", [False, True], ids=["tau8", "exact_max"])
def test_pair64_row_max_rising_across_tiles(exact):
    """Keys scaled up along the sequence, so each row's max rises tile after
    tile; in exact-max mode O is rescaled on most tiles."""
    q, k, v = inputs.make_qkv(1, 4, 1100, 1100, 128, "fp16", 35, qk_mult=2.0)
    ramp = 1.0 + 3.0 * torch.arange(k.shape[2], dtype=torch.float32) / k.shape[2]
    k = (k.float() * ramp[None, None, :, None]).to(k.dtype)
    f = P64 | (fa.FA_FLAG_EXACT_MAX if exact else 0)
    o, lse = run_kernel(q, k, v, False, flags=f)
    _assert(check(q, k, v, o, lse, False, "fp16"))
    o2, l2 = run_kernel(q, k, v, False, flags=f | fa.FA_FLAG_ALWAYS_RESCALE)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_pair64_watchdog_reports_timeout_and_context_survives():
    q, k, v = inputs.make_qkv(1, 2, 512, 512, 128, "bf16", 36)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)
    try:
        fa.fa_fwd_ex(dq, dk, dv, flags=P64 | fa.FA_FLAG_TEST_STALL)
        assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_device_status() == fa.FA_OK
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = run_kernel(q, k, v, False, flags=P64)
    _assert(check(q, k, v, o, lse, False, "bf16"))
