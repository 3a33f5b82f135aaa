"""Parity of the three-stage D = 64 prefill kernel (FA_FLAG_D64_THREE_STAGE:
384-row items of three 128-row stages, 96-key tiles) with the fp64 oracle,
through the C ABI.  Gate: oracle/gate.py."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_and_check, run_kernel, sample_rows

pytestmark = pytest.mark.gpu

X3 = fa.FA_FLAG_D64_THREE_STAGE


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _assert(r):
    assert r.passed, str(r)


CASES = [  # B, H, Sq, Skv, dtype, causal
    (1, 1, 2, 2, "bf16", True),        # one item, almost all rows padding
    (1, 1, 96, 96, "fp16", False),     # one key tile exactly
    (1, 1, 97, 97, "bf16", True),      # a ragged second tile
    (1, 2, 129, 129, "bf16", True),    # stage 2 past Sq, stage 1 one row
    (1, 1, 256, 300, "fp16", False),   # stage 2 past Sq
    (1, 1, 383, 383, "bf16", True),
    (1, 1, 384, 384, "bf16", False),   # one full item
    (1, 1, 385, 385, "fp16", True),    # two items, the second one row
    (2, 3, 1000, 1000, "bf16", True),
    (1, 1, 100, 300, "fp16", True),    # Sq < Skv (bottom-right diagonal)
    (1, 1, 300, 100, "bf16", True),    # Sq > Skv: rows without a visible key
    (1, 1, 600, 40, "bf16", False),    # fewer keys than one tile
    (1, 1, 800, 129, "fp16", True),
    (2, 8, 1024, 1024, "bf16", False),
    (2, 8, 1024, 1024, "bf16", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_d64x3_edge_shapes(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 64, dt, causal, 41, qk_mult=2.0, flags=X3))


# more items than SMs: every CTA takes several items in turn
PERSISTENT = [
    (4, 48, 600, 129, "bf16", True),
    (8, 32, 300, 300, "bf16", False),
    (1, 64, 1024, 128, "fp16", True),
    (4, 16, 2048, 2048, "bf16", True),
    (2, 16, 2048, 2048, "fp16", False),
]


@pytest.mark.parametrize("case", PERSISTENT, ids=lambda c: "x".join(map(str, c)))
def test_d64x3_persistent_item_sequences(case):
    B, H, Sq, Skv, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, 64, dt, causal, 42, flags=X3))


@pytest.mark.parametrize("name", ["sweep_S4096_D64_bf16_full", "sweep_S4096_D64_bf16_causal",
                                  "sweep_S16384_D64_fp16_causal"])
def test_d64x3_sweep_sampled_rows(name):
    w = inputs.BY_NAME[name]
    rows = sample_rows(w.B, w.H, w.Sq, per_head=24, extra=256, seed=9)
    assert rows.size >= 512
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed,
                          rows=rows, flags=X3))


def test_d64x3_repeat_and_switches_bitwise_identical():
    """Repeats, the plain item order and rescaling on every tile give the
    same bits."""
    q, k, v = inputs.make_qkv(4, 16, 1500, 1500, 64, "bf16", 43, 4.0)
    o1, l1 = run_kernel(q, k, v, True, flags=X3)
    o2, l2 = run_kernel(q, k, v, True, flags=X3)
    o3, l3 = run_kernel(q, k, v, True, flags=X3 | fa.FA_FLAG_NO_LPT)
    o4, l4 = run_kernel(q, k, v, True, flags=X3 | fa.FA_FLAG_ALWAYS_RESCALE)
    for o, l in ((o2, l2), (o3, l3), (o4, l4)):
        assert torch.equal(o, o1) and torch.equal(l, l1)


@pytest.mark.parametrize("scale", [1.0, 1e-3], ids=["sharp", "flat"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_d64x3_extreme_scales(scale, causal):
    q, k, v = inputs.make_qkv(1, 4, 1500, 1500, 64, "bf16", 44)
    v = v * 0.25
    o, lse = run_kernel(q, k, v, causal, flags=X3, scale=scale)
    _assert(check(q, k, v, o, lse, causal, "bf16", scale=scale))


@pytest.mark.parametrize("exact", [False, True], ids=["tau8", "exact_max"])
def test_d64x3_row_max_rising_across_tiles(exact):
    q, k, v = inputs.make_qkv(1, 4, 1100, 1100, 64, "fp16", 45, qk_mult=2.0)
    ramp = 1.0 + 3.0 * torch.arange(k.shape[2], dtype=torch.float32) / k.shape[2]
    k = (k.float() * ramp[None, None, :, None]).to(k.dtype)
    f = X3 | (fa.FA_FLAG_EXACT_MAX if exact else 0)
    o, lse = run_kernel(q, k, v, False, flags=f)
    _assert(check(q, k, v, o, lse, False, "fp16"))
    o2, l2 = run_kernel(q, k, v, False, flags=f | fa.FA_FLAG_ALWAYS_RESCALE)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_d64x3_overlapped_calls_match_plain_calls():
    q, k, v = (t.cuda() for t in inputs.make_qkv(4, 16, 2048, 2048, 64, "bf16", 46))
    ref_o, ref_l = fa.fa_fwd_ex(q, k, v, causal=True, flags=X3)
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    for _ in range(20):
        fa.fa_fwd_ex(q, k, v, causal=True, flags=X3 | fa.FA_FLAG_OVERLAP_PREVIOUS, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_d64x3_flag_ignored_where_it_does_not_apply():
    """D = 128 and an explicit key split run the other kernels."""
    _assert(run_and_check(1, 2, 300, 300, 128, "bf16", True, 47, flags=X3))
    q, k, v = inputs.make_qkv(1, 2, 256, 2048, 64, "bf16", 48)
    need = fa.fa_workspace_bytes(1, 2, 256, 2048, 64, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = run_kernel(q, k, v, True, flags=X3, num_splits=4, workspace=ws)
    _assert(check(q, k, v, o, lse, True, "bf16"))


def test_d64x3_watchdog_reports_timeout_and_context_survives():
    q, k, v = inputs.make_qkv(1, 2, 512, 512, 64, "bf16", 49)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)
    try:
        fa.fa_fwd_ex(dq, dk, dv, flags=X3 | fa.FA_FLAG_TEST_STALL)
        assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_device_status() == fa.FA_OK
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = run_kernel(q, k, v, False, flags=X3)
    _assert(check(q, k, v, o, lse, False, "bf16"))
